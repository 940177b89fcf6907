"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (bulk tq_quantize_kv of the whole context, then
tq_decode_attention over every sequence and head with one workspace).

The oracle cannot redo a whole full-size call in seconds, so it recomputes
sampled (sequence, kv-head) pairs one by one from the same seeded inputs:
their packed codes (bit-exact but for the boundary band) and the attention
output of the kv-head's query heads (2e-3 relative L2).
"""

import numpy as np
import pytest

import oracle as O
from gpu_helpers import binding, rel_l2_per_head, to64

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def B():
    return binding()


def _layer_cache(B, w, cfg, tables, layer, seq, device):
    """Seeded K/V of one layer on the GPU, bulk-quantized into planes, plus the
    bf16 window ring of every sequence."""
    import torch
    from kv_cache_quantization_random_gb300 import workloads as WL
    K, V = WL.make_kv(w, layer=layer, device=device)
    Wn = w.window
    Tmax = int(seq.max())
    nq = max(Tmax - Wn, 0)
    kp = B.Planes(cfg, layer, 0, w.batch, w.n_kv_heads, max(nq, 1), device)
    vp = B.Planes(cfg, layer, 1, w.batch, w.n_kv_heads, max(nq, 1), device)
    if nq:
        B.tq_quantize_kv(cfg, tables, layer, 0, K[:, :, :nq], kp)
        B.tq_quantize_kv(cfg, tables, layer, 1, V[:, :, :nq], vp)
    kw = vw = None
    if Wn:
        kw = torch.zeros(w.batch, w.n_kv_heads, Wn, w.head_dim, dtype=torch.bfloat16, device=device)
        vw = torch.zeros_like(kw)
        for b in range(w.batch):
            T = int(seq[b])
            t = torch.arange(max(T - Wn, 0), T, device=device)
            kw[b, :, t % Wn] = K[b, :, t]
            vw[b, :, t % Wn] = V[b, :, t]
    return K, V, kp, vp, kw, vw


def _check_samples(B, w, cfg, layer, K, V, kp, vp, q, out, seq, samples):
    """Oracle quantize + decode of each sampled (b, kv-head) against the GPU."""
    kb, vb, mode = B.tq_layer_spec_get(cfg, layer)
    seed = w.codec_seed
    ck, bk = O.codebook_fp32(kb, w.head_dim)
    cv, bv = O.codebook_fp32(vb, w.head_dim)
    sk = O.rotation_signs(seed, layer, 0, w.head_dim)
    sv = O.rotation_signs(seed, layer, 1, w.head_dim)
    g = w.group
    Wn = w.window
    worst = 0.0
    for b, h in samples:
        T = int(seq[b])
        nq = max(T - Wn, 0)
        K64 = to64(K[b:b + 1, h:h + 1, :T])
        V64 = to64(V[b:b + 1, h:h + 1, :T])
        qk = O.quantize_vectors(K64[:, :, :nq], ck, bk, sk)
        qv = O.quantize_vectors(V64[:, :, :nq], cv, bv, sv)
        # codes: every row up to 65,536 rows, else an evenly strided subset
        rows = np.arange(nq)[::max(1, nq // 65536)]
        for planes, oq, bits, b32 in ((kp, qk, kb, bk), (vp, qv, vb, bv)):
            gpu = O.unpack_codes(planes.codes_view()[b, h].cpu().numpy()[rows], bits, w.head_dim)
            ref_codes = oq["codes"][0, 0][rows]
            diff = gpu != ref_codes
            if diff.any():
                band = O.near_boundary(oq["y"][0, 0][rows][diff], b32, w.head_dim)
                assert band.all(), int((~band).sum())
                assert np.abs(gpu[diff] - ref_codes[diff]).max() <= 1
        qjl = None
        if mode == B.TQ_MODE_MSE_QJL:
            S = O.qjl_matrix(seed, layer, w.qjl_m, w.head_dim)
            r = O.qjl_residual(qk["y"], qk["codes"], qk["norm64"], ck)
            bits, gamma, _ = O.qjl_sketch(r, S)
            qjl = dict(bits=bits, gamma=gamma, S=S)
        kw = vw = None
        if Wn:
            kw = np.zeros((1, 1, Wn, w.head_dim))
            vw = np.zeros_like(kw)
            for t in range(nq, T):
                kw[0, 0, t % Wn] = K64[0, 0, t]
                vw[0, 0, t % Wn] = V64[0, 0, t]
        qs = to64(q[b:b + 1, h * g:(h + 1) * g])
        ref = O.decode_attention(qs, qk["codes"], qk["norms"], qv["codes"], qv["norms"], ck, cv,
                                 sk, sv, [T], w.softmax_scale, window=Wn, k_win=kw, v_win=vw,
                                 qjl=qjl)
        got = to64(out[b:b + 1, h * g:(h + 1) * g])
        rel = rel_l2_per_head(got, ref).max()
        worst = max(worst, float(rel))
        assert rel < TOL, (b, h, rel)
    return worst


def _decode(B, w, cfg, tables, layer, kp, vp, kw, vw, seq, device):
    import torch
    from kv_cache_quantization_random_gb300 import workloads as WL
    q = WL.make_q(w, layer=layer, device=device)
    Tmax = int(seq.max())
    out = torch.full((w.batch, w.n_q_heads, w.head_dim), float("nan"), device=device)
    ws = B.new_workspace(cfg, w.batch, w.n_q_heads, w.n_kv_heads, Tmax, device)
    seq_t = torch.tensor(seq, dtype=torch.int32, device=device)
    B.tq_decode_attention(cfg, tables, layer, q, w.softmax_scale, kp, vp, seq_t, Tmax, out, ws,
                          k_win=kw, v_win=vw)
    torch.cuda.synchronize()
    assert B.tq_get_device_error() == B.TQ_OK
    assert torch.isfinite(out).all()
    return q, out


@pytest.mark.parametrize("name", ["llama8b_32k", "qjl_b16_8k", "long_1m"])
def test_full_size_quantize_and_decode(B, name):
    import torch
    from kv_cache_quantization_random_gb300 import workloads as WL
    w = WL.get(name)
    dev = torch.device("cuda", 0)
    cfg = B.Config(k_bits=w.k_bits, v_bits=w.v_bits, residual_window=w.window, seed=w.codec_seed,
                   k_mode=B.TQ_MODE_MSE_QJL if w.k_qjl else B.TQ_MODE_MSE, qjl_m=w.qjl_m)
    tables = B.device_tables(cfg, dev)
    seq = WL.seq_lens(w)
    K, V, kp, vp, kw, vw = _layer_cache(B, w, cfg, tables, 0, seq, dev)
    q, out = _decode(B, w, cfg, tables, 0, kp, vp, kw, vw, seq, dev)
    samples = [(0, 0), (w.batch - 1, w.n_kv_heads - 1)]
    if name == "long_1m":
        samples = [(0, 3)]              # one kv-head of the 1M-token sequence
    _check_samples(B, w, cfg, 0, K, V, kp, vp, q, out, seq, samples)


def test_serving_36_layers_full_batch(B):
    """The 36-layer serving stack at full batch (64 ragged sequences of 4K-16K
    tokens): protected 8-bit layers and K4/V2 layers, sampled per layer."""
    import torch
    from kv_cache_quantization_random_gb300 import workloads as WL
    w = WL.get("serving_36l")
    dev = torch.device("cuda", 0)
    cfg = B.Config(n_layers=w.n_layers, k_bits=w.k_bits, v_bits=w.v_bits,
                   n_protect_first=w.protect_first, n_protect_last=w.protect_last,
                   residual_window=w.window, seed=w.codec_seed)
    tables = B.device_tables(cfg, dev)
    seq = WL.seq_lens(w)
    shortest, longest = int(np.argmin(seq)), int(np.argmax(seq))
    for layer in (0, 4, 35):
        K, V, kp, vp, kw, vw = _layer_cache(B, w, cfg, tables, layer, seq, dev)
        q, out = _decode(B, w, cfg, tables, layer, kp, vp, kw, vw, seq, dev)
        samples = [(shortest, 0), (longest, w.n_kv_heads - 1), (w.batch // 2, 3)]
        _check_samples(B, w, cfg, layer, K, V, kp, vp, q, out, seq, samples)
        del K, V, kp, vp
        torch.cuda.empty_cache()
