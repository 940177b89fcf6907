"""The allocation-free decode entry point (tq_decode_attention_noalloc).

Some callers cannot hand the library a workspace: a plugin inside a serving
engine that owns every device allocation and passes only tensor pointers, or
a latency-bound decode loop that must not call the CUDA allocator (cudaMalloc
can synchronize the whole device).  This entry point keeps the decode scratch
in a fixed device array inside the library instead.

The GPU test runs two calls in a row with different shapes (so what the first
call leaves in the shared array must not leak into the second).  Each output
must be bit-identical to tq_decode_attention with a caller workspace (the same
kernel runs the same split plan) and within the decode tolerance of the oracle,
run on the oracle's own quantization of the same seeded inputs.  A host test
checks that an oversized problem is refused before anything is launched.  The
file is named so that pytest collects it last.
"""

import ctypes as C

import numpy as np
import pytest

from gpu_helpers import rel_l2_per_head

TOL = 2e-3


@pytest.mark.gpu
def test_noalloc_decode_matches_workspace_decode_and_oracle_on_two_calls():
    import torch
    from gpu_helpers import binding
    from test_gpu_decode import _decode_case
    B = binding()
    cases = [
        dict(batch=2, hq=8, hkv=2, seq=[1500, 333], kb=4, vb=2, W=16, data_seed=21),
        dict(batch=3, hq=16, hkv=2, seq=[17, 900, 500], kb=3, vb=3, W=32, data_seed=22),
    ]
    for case in cases:      # two calls in a row, different shapes
        ws_out, ref, c = _decode_case(B, **case)
        got = torch.full((case["batch"], case["hq"], 128), float("nan"), device="cuda")
        B.tq_decode_attention_noalloc(c["cfg"], c["tables"], 0, c["q"].cuda(), c["scale"],
                                      c["kp"], c["vp"], c["seq_t"], c["Tmax"], got,
                                      k_win=c["kw"], v_win=c["vw"])
        torch.cuda.synchronize()
        assert B.tq_get_device_error() == B.TQ_OK
        g = got.double().cpu().numpy()
        assert np.array_equal(g, ws_out)
        assert rel_l2_per_head(g, ref).max() < TOL


def test_noalloc_rejects_problems_larger_than_its_array():
    """Host-side size check: the call must refuse before any memset or launch,
    so it never touches the (tiny) buffers it is given."""
    from conftest import has_gpu
    from kv_cache_quantization_random_gb300 import binding as B
    from kv_cache_quantization_random_gb300 import build
    if not has_gpu():
        build.build()
    lib = B.load(build_if_missing=True)
    cfg = B.Config(residual_window=128)
    batch, hq, hkv, T = 256, 64, 8, 1 << 20
    assert B.tq_workspace_bytes(cfg, batch, hq, hkv, T) > B.NOALLOC_MAX_BYTES
    if has_gpu():
        import torch
        buf = torch.zeros(64, dtype=torch.float32, device="cuda")     # 256 bytes, never read
        p = buf.data_ptr()
    else:
        p = 4096                                                       # placeholder, never read
    planes = B.tq_planes(p, p, None, None, T)
    rc = lib.tq_decode_attention_noalloc(C.byref(cfg.c()), p, 0, p, 0, 1.0, batch, hq, hkv,
                                         planes, planes, p, p, p, T, p, None)
    assert rc == B.TQ_ERR_BUFFER_TOO_SMALL
