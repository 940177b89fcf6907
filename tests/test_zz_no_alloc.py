"""The allocation-free decode entry point (tq_decode_attention_noalloc).

Callers such as a plugin inside a serving engine that owns all device memory,
or a latency-bound decode loop that must not call the CUDA allocator, cannot
pass a workspace; this entry point keeps the decode scratch in a fixed device
array inside the library instead.  These tests check that it gives the same
attention output as tq_decode_attention with a caller workspace, on two calls
in a row with different problem sizes (so leftovers of the first call in the
shared array must not leak into the second), and that an oversized problem is
rejected before anything runs.  The file is named so that pytest collects it
last.
"""

import ctypes as C

import numpy as np
import pytest

TOL = 2e-3


def _rel_l2(a, b):
    num = np.linalg.norm(a - b, axis=-1)
    den = np.linalg.norm(b, axis=-1)
    return np.where(den > 0, num / np.maximum(den, 1e-300), num)


def _cache(B, torch, batch, hq, hkv, T, W, seed):
    from kv_cache_quantization_random_gb300 import workloads as WL
    w = WL.scaled(WL.get("llama8b_32k"), batch=batch, n_q_heads=hq, n_kv_heads=hkv, context=T,
                  window=W, data_seed=seed)
    K, V = WL.make_kv(w)
    nq = T - W
    cfg = B.Config(k_bits=4, v_bits=2, residual_window=W, seed=seed)
    tables = B.device_tables(cfg)
    kp = B.Planes(cfg, 0, 0, batch, hkv, nq)
    vp = B.Planes(cfg, 0, 1, batch, hkv, nq)
    B.tq_quantize_kv(cfg, tables, 0, 0, K[:, :, :nq].cuda(), kp)
    B.tq_quantize_kv(cfg, tables, 0, 1, V[:, :, :nq].cuda(), vp)
    kw = torch.empty(batch, hkv, W, 128, dtype=torch.bfloat16)
    vw = torch.empty_like(kw)
    for t in range(nq, T):
        kw[:, :, t % W] = K[:, :, t]
        vw[:, :, t % W] = V[:, :, t]
    return dict(w=w, cfg=cfg, tables=tables, kp=kp, vp=vp, kw=kw.cuda(), vw=vw.cuda(),
                q=WL.make_q(w).cuda())


@pytest.mark.gpu
def test_noalloc_decode_matches_workspace_decode_on_two_calls():
    import torch
    from kv_cache_quantization_random_gb300 import binding as B
    B.load(build_if_missing=True)
    cases = [
        dict(batch=2, hq=8, hkv=2, T=1500, W=16, seed=21, seq=[1500, 333]),
        dict(batch=3, hq=16, hkv=2, T=900, W=32, seed=22, seq=[17, 900, 500]),
    ]
    for case in cases:      # two calls in a row, different shapes
        c = _cache(B, torch, case["batch"], case["hq"], case["hkv"], case["T"], case["W"],
                   case["seed"])
        seq = torch.tensor(case["seq"], dtype=torch.int32, device="cuda")
        Tmax = max(case["seq"])
        ref = torch.empty(case["batch"], case["hq"], 128, device="cuda")
        ws = B.new_workspace(c["cfg"], case["batch"], case["hq"], case["hkv"], Tmax)
        B.tq_decode_attention(c["cfg"], c["tables"], 0, c["q"], c["w"].softmax_scale, c["kp"],
                              c["vp"], seq, Tmax, ref, ws, k_win=c["kw"], v_win=c["vw"])
        got = torch.full_like(ref, float("nan"))
        B.tq_decode_attention_noalloc(c["cfg"], c["tables"], 0, c["q"], c["w"].softmax_scale,
                                      c["kp"], c["vp"], seq, Tmax, got, k_win=c["kw"],
                                      v_win=c["vw"])
        torch.cuda.synchronize()
        assert B.tq_get_device_error() == B.TQ_OK
        r = ref.double().cpu().numpy()
        g = got.double().cpu().numpy()
        assert np.all(np.isfinite(g))
        assert _rel_l2(g, r).max() < TOL


def test_noalloc_rejects_problems_larger_than_its_array():
    """Host-side size check (runs without a GPU: it must refuse before any launch)."""
    from conftest import has_gpu
    if has_gpu():
        pytest.skip("uses placeholder pointers, which only a machine without a GPU may see")
    from kv_cache_quantization_random_gb300 import binding as B
    from kv_cache_quantization_random_gb300 import build
    build.build()
    lib = B.load()
    cfg = B.Config(residual_window=128)
    batch, hq, hkv, T = 256, 64, 8, 1 << 20
    assert B.tq_workspace_bytes(cfg, batch, hq, hkv, T) > B.NOALLOC_MAX_BYTES
    planes = B.tq_planes(4096, 8192, None, None, T)
    rc = lib.tq_decode_attention_noalloc(C.byref(cfg.c()), 4096, 0, 16384, 0, 1.0, batch, hq,
                                         hkv, planes, planes, 32768, 32768, 20480, T, 65536, None)
    assert rc == 7          # TQ_ERR_BUFFER_TOO_SMALL
