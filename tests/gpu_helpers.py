"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same seeded inputs, compare."""

import math

import numpy as np

import oracle as O


def binding():
    from kv_cache_quantization_random_gb300 import binding as B
    B.load(build_if_missing=True)
    return B


def to64(t):
    """Exact fp64 copy of a torch tensor (bf16 / fp32)."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def oracle_codec(bits, d=128):
    return O.codebook_fp32(bits, d)


def oracle_codebook(bits, d=128, density=0):
    """fp32 codebook of the oracle: N(0, 1/d) (density 0) or sphere (1)."""
    return O.codebook_sphere_fp32(bits, d) if density == 1 else O.codebook_fp32(bits, d)


def oracle_quantize(X64, bits, seed, layer, kind, d=128, density=0):
    c32, b32 = oracle_codebook(bits, d, density)
    s = O.rotation_signs(seed, layer, kind, d)
    q = O.quantize_vectors(X64, c32, b32, s)
    q["packed"] = O.pack_codes(q["codes"], bits)
    q["c32"], q["b32"], q["signs"] = c32, b32, s
    return q


def compare_codes(gpu_packed, oq, bits, d=128):
    """Packed codes must be bit-exact, except coordinates within 1e-6 relative
    of a decision boundary, which may differ by one code.  Returns the number of
    such coordinates."""
    gpu_codes = O.unpack_codes(gpu_packed, bits, d)
    diff = gpu_codes != oq["codes"]
    if diff.any():
        band = O.near_boundary(oq["y"], oq["b32"], d, rel=1e-6)
        bad = diff & ~band
        assert not bad.any(), f"{int(bad.sum())} code mismatches outside the boundary band"
        assert np.abs(gpu_codes - oq["codes"])[diff].max() <= 1
    else:
        assert np.array_equal(gpu_packed, oq["packed"])
    return int(diff.sum())


def compare_norms(gpu, oracle32, rel=1e-6):
    g = np.asarray(gpu, dtype=np.float64)
    o = np.asarray(oracle32, dtype=np.float64)
    err = np.abs(g - o)
    assert np.all(err <= rel * np.abs(o) + 1e-30), float((err / np.maximum(np.abs(o), 1e-30)).max())


def rel_l2_per_head(out, ref):
    num = np.linalg.norm(out - ref, axis=-1)
    den = np.linalg.norm(ref, axis=-1)
    return np.where(den > 0, num / np.maximum(den, 1e-300), num)


def upload_oracle_planes(B, planes, oq, layer_rows=None):
    """Write the oracle's packed codes / fp32 norms into GPU planes
    (rows [0, T) of every (sequence, head))."""
    import torch
    Bsz, H, T = oq["codes"].shape[:3]
    cv = planes.codes_view()
    cv[:, :, :T].copy_(torch.from_numpy(np.ascontiguousarray(oq["packed"])))
    planes.norms_view()[:, :, :T].copy_(torch.from_numpy(np.ascontiguousarray(oq["norms"])))


def oracle_qjl(oq, seed, layer, m=128, d=128):
    S = O.qjl_matrix(seed, layer, m, d)
    r = O.qjl_residual(oq["y"], oq["codes"], oq["norm64"], oq["c32"])
    bits, gamma, z = O.qjl_sketch(r, S)
    return dict(S=S, bits=bits, gamma=gamma, z=z, packed=O.pack_bits(bits), r=r)


def oq_slice(oq, idx):
    """The oracle result restricted to an index expression over its leading axes."""
    return dict(codes=oq["codes"][idx], y=oq["y"][idx], packed=oq["packed"][idx],
                norms=oq["norms"][idx], b32=oq["b32"], c32=oq["c32"], signs=oq["signs"])
