"""Seeded synthetic workloads: shapes, sizes and value distributions only.

This module holds none of the codec's arithmetic.  It is the one module that
both the CUDA path's tests and benchmark and the CPU oracle's inputs come from.

The five workloads mirror the shapes on the TurboQuant pages:

* ``single_head_1k``  one head, d = 128, 1024 tokens, fp32 K/V ~ N(0,1) with 4
  outlier channels x20, 3-bit keys and values, query N(0,1)/sqrt(d) (already
  scaled, so the softmax scale is 1).
* ``llama8b_32k``  Llama-3-8B-shaped decode layer: batch 1, 32 query / 8 KV
  heads, 32768 tokens, bf16; keys with log-normal(0,1) per-channel sigma, 6
  outlier channels (5 % of 128) x20, rescaled to a mean key norm of about 170;
  values N(0, 0.25^2) (norm about 3); K4/V2, residual window of 128 tokens.
  The key/value norm gap is the one the write-up measured on Qwen2.5 caches
  ("윈도우용 터보퀀트(TurboQuant) 구현을 개선하다", finding 2).
* ``qjl_b16_8k``  batch 16, 32/8 heads, 8192 tokens, keys 2-bit + 1-bit QJL
  sketch (m = 128), values 3-bit, no window.
* ``sign_b16_8k``  the same shapes and inputs with the keys' 1-bit residual
  term stored as Direct Sign (128 residual signs + scale) instead of QJL.
* ``long_1m``  batch 1, 64/8 heads, 1,048,576 tokens, K3/V3, window 256,
  streaming quantize in 4096-token chunks.
* ``serving_36l``  36 layers, layers 0-3 and 32-35 at 8 bits, the rest K4/V2;
  batch 64, 32/8 heads, contexts uniform in [4096, 16384], 64 new tokens per
  sequence per step.
The QJL, Direct Sign, long-context and serving workloads draw their keys and
values from the first workload's distributions (N(0,1) with 4 outlier channels
x20, keys and values alike), in bf16, with a query N(0,1) and softmax scale
1/sqrt(d).  ``with_llama_kv`` gives the same shapes with the Llama-shaped
key/value distributions instead (a bench option).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional, Tuple

import numpy as np

__all__ = ["Workload", "WORKLOADS", "get", "seq_lens", "kv_params", "make_kv", "make_q",
           "scaled", "with_llama_kv"]


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    context: int                       # tokens per sequence (max when ragged)
    k_bits: int
    v_bits: int
    k_qjl: bool = False
    k_sign: bool = False               # keys with the Direct Sign residual
    qjl_m: int = 128
    window: int = 0
    n_layers: int = 1
    protect_first: int = 0
    protect_last: int = 0
    protect_bits: int = 8
    in_dtype: str = "bf16"             # "bf16" | "fp32"
    dist: str = "llama"                # "gauss_outlier" | "llama"
    n_outliers: int = 6
    outlier_gain: float = 20.0
    key_norm: float = 170.0
    value_sigma: float = 0.25
    query_prescaled: bool = False      # q ~ N(0,1)/sqrt(d) and softmax scale 1
    ragged: Optional[Tuple[int, int]] = None
    new_tokens: int = 1                # tokens appended per decode step
    data_seed: int = 1000
    codec_seed: int = 0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def softmax_scale(self) -> float:
        return 1.0 if self.query_prescaled else 1.0 / math.sqrt(self.head_dim)


WORKLOADS = {
    "single_head_1k": Workload(
        name="single_head_1k", batch=1, n_q_heads=1, n_kv_heads=1, head_dim=128,
        context=1024, k_bits=3, v_bits=3, in_dtype="fp32", dist="gauss_outlier",
        n_outliers=4, query_prescaled=True, data_seed=1000),
    "llama8b_32k": Workload(
        name="llama8b_32k", batch=1, n_q_heads=32, n_kv_heads=8, head_dim=128,
        context=32768, k_bits=4, v_bits=2, window=128, data_seed=1001),
    "qjl_b16_8k": Workload(
        name="qjl_b16_8k", batch=16, n_q_heads=32, n_kv_heads=8, head_dim=128,
        context=8192, k_bits=2, v_bits=3, k_qjl=True, qjl_m=128, data_seed=1002,
        dist="gauss_outlier", n_outliers=4),
    "sign_b16_8k": Workload(
        name="sign_b16_8k", batch=16, n_q_heads=32, n_kv_heads=8, head_dim=128,
        context=8192, k_bits=2, v_bits=3, k_sign=True, data_seed=1002,
        dist="gauss_outlier", n_outliers=4),
    "long_1m": Workload(
        name="long_1m", batch=1, n_q_heads=64, n_kv_heads=8, head_dim=128,
        context=1048576, k_bits=3, v_bits=3, window=256, new_tokens=4096,
        data_seed=1003,
        dist="gauss_outlier", n_outliers=4),
    "serving_36l": Workload(
        name="serving_36l", batch=64, n_q_heads=32, n_kv_heads=8, head_dim=128,
        context=16384, k_bits=4, v_bits=2, n_layers=36, protect_first=4,
        protect_last=4, ragged=(4096, 16384), new_tokens=64, data_seed=1004,
        dist="gauss_outlier", n_outliers=4),
}


def get(name: str) -> Workload:
    return WORKLOADS[name]


def with_llama_kv(w: Workload) -> Workload:
    """The same shapes with the Llama-shaped key/value distributions
    (log-normal key channels, 6 outliers, mean key norm 170, values
    N(0, 0.25^2))."""
    return replace(w, dist="llama", n_outliers=6)


def scaled(w: Workload, **kw) -> Workload:
    """The same workload with some sizes changed (small parity cases)."""
    return replace(w, **kw)


def seq_lens(w: Workload) -> np.ndarray:
    """Tokens per sequence (window included), int32 [batch]."""
    if w.ragged is None:
        return np.full(w.batch, w.context, dtype=np.int32)
    rng = np.random.default_rng(w.data_seed + 17)
    lo, hi = w.ragged
    return rng.integers(lo, hi + 1, size=w.batch).astype(np.int32)


def kv_params(w: Workload, layer: int = 0):
    """Per-(kv-head, channel) key scale and value scale, [Hkv, d] float64.

    llama: sigma_c = exp(N(0,1)); n_outliers channels (without replacement)
    x outlier_gain; the head is then rescaled so that the mean key norm is
    key_norm.  gauss_outlier: unit sigma with outliers, applied to
    keys and values alike.
    """
    rng = np.random.default_rng([w.data_seed, layer, 7])
    H, d = w.n_kv_heads, w.head_dim
    ks = np.empty((H, d))
    vs = np.empty((H, d))
    for h in range(H):
        out = rng.choice(d, size=w.n_outliers, replace=False)
        if w.dist == "llama":
            sig = np.exp(rng.standard_normal(d))
            sig[out] *= w.outlier_gain
            # rescale so that the mean key norm is key_norm: the norm of
            # sigma * z has no closed-form mean, so measure it on a fixed
            # seeded sample of 4096 vectors
            probe = np.random.default_rng([w.data_seed, layer, h, 11]).standard_normal((4096, d))
            sig *= w.key_norm / np.mean(np.linalg.norm(probe * sig, axis=1))
            ks[h] = sig
            vs[h] = w.value_sigma
        elif w.dist == "gauss_outlier":
            sig = np.ones(d)
            sig[out] *= w.outlier_gain
            ks[h] = sig
            vs[h] = sig
        else:
            raise ValueError(w.dist)
    return ks, vs


def _torch_dtype(w: Workload):
    import torch
    return torch.float32 if w.in_dtype == "fp32" else torch.bfloat16


def make_kv(w: Workload, layer: int = 0, device="cpu", tokens: Optional[int] = None,
            batch: Optional[int] = None, token_offset: int = 0):
    """K and V as torch tensors [B, Hkv, T, d] in the workload's input dtype.

    The noise comes from a torch generator seeded by (data_seed, layer,
    token_offset), on ``device``; drawing the same slice twice on the same
    device gives the same tensors.
    """
    import torch
    T = w.context if tokens is None else tokens
    B = w.batch if batch is None else batch
    ks, vs = kv_params(w, layer)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(w.data_seed) * 1_000_003 + layer * 7919 + token_offset)
    shape = (B, w.n_kv_heads, T, w.head_dim)
    K = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    K.mul_(torch.as_tensor(ks, dtype=torch.float32, device=device)[None, :, None, :])
    V = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    V.mul_(torch.as_tensor(vs, dtype=torch.float32, device=device)[None, :, None, :])
    dt = _torch_dtype(w)
    return K.to(dt), V.to(dt)


def make_q(w: Workload, layer: int = 0, device="cpu", step: int = 0):
    """Decode queries [B, Hq, d]: N(0,1), or N(0,1)/sqrt(d) when prescaled."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(w.data_seed) * 999_983 + layer * 31 + step)
    q = torch.randn((w.batch, w.n_q_heads, w.head_dim), generator=gen, device=device,
                    dtype=torch.float32)
    if w.query_prescaled:
        q.mul_(1.0 / math.sqrt(w.head_dim))
    return q.to(_torch_dtype(w))
