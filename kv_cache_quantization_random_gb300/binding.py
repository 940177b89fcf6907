"""Thin Python binding of the TurboQuant C ABI (include/tq.h).

Argument marshalling only: every step of the path runs in the CUDA library.
PyTorch provides device memory and streams.  The functions carry the C names
(``tq_quantize_kv`` ...) and take torch tensors where the C call takes device
pointers.  There is no CPU fallback: if ``libtq.so`` is missing, loading fails
with an error that says how to build it.
"""

from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

from . import build as _build

TQ_OK = 0
TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_ALIGNMENT, TQ_ERR_CUDA = 1, 2, 3, 4
TQ_ERR_DEVICE_TIMEOUT, TQ_ERR_DEVICE_BOUNDS, TQ_ERR_BUFFER_TOO_SMALL = 5, 6, 7
TQ_ERR_NAMES = {
    0: "TQ_OK", 1: "TQ_ERR_INVALID_ARG", 2: "TQ_ERR_UNSUPPORTED", 3: "TQ_ERR_ALIGNMENT",
    4: "TQ_ERR_CUDA", 5: "TQ_ERR_DEVICE_TIMEOUT", 6: "TQ_ERR_DEVICE_BOUNDS",
    7: "TQ_ERR_BUFFER_TOO_SMALL",
}
TQ_MODE_MSE, TQ_MODE_MSE_QJL, TQ_MODE_MSE_SIGN = 0, 1, 2
TQ_DENSITY_GAUSSIAN, TQ_DENSITY_SPHERE_BETA = 0, 1
TQ_BF16, TQ_F32 = 0, 1
TQ_KIND_K, TQ_KIND_V = 0, 1

# every symbol include/tq.h declares
EXPORTED = [
    "tq_version", "tq_status_string", "tq_layer_spec_get", "tq_make_codebook", "tq_make_signs",
    "tq_make_qjl_matrix", "tq_tables_bytes", "tq_build_tables", "tq_plane_bytes",
    "tq_workspace_bytes", "tq_workspace_init", "tq_quantize_kv", "tq_append_kv",
    "tq_dequantize", "tq_decode_attention", "tq_get_device_error", "tq_set_wait_limit",
    "tq_set_fault_injection", "tq_decode_attention_noalloc", "tq_decode_attention_multi",
    "tq_decode_step", "tq_decode_step_launches",
]


class TQError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {TQ_ERR_NAMES.get(status, status)}")
        self.status = status


class tq_config(C.Structure):
    _fields_ = [("head_dim", C.c_int32), ("n_layers", C.c_int32), ("k_bits", C.c_int32),
                ("v_bits", C.c_int32), ("k_mode", C.c_int32), ("qjl_m", C.c_int32),
                ("n_protect_first", C.c_int32), ("n_protect_last", C.c_int32),
                ("protect_bits", C.c_int32), ("residual_window", C.c_int32),
                ("density", C.c_int32), ("sparse_v", C.c_int32), ("seed", C.c_uint64)]


class tq_layer_spec(C.Structure):
    _fields_ = [("k_bits", C.c_int32), ("v_bits", C.c_int32), ("k_mode", C.c_int32)]


class tq_planes(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("norms", C.c_void_p), ("qjl_signs", C.c_void_p),
                ("qjl_rnorm", C.c_void_p), ("capacity", C.c_int64)]


_LIB = None


def lib_path() -> str:
    """The library this process loads: libtq.so, or with TQ_LIB_VARIANT=debug
    the bounds-checked libtq_debug.so."""
    return _build.lib_path()


def load(build_if_missing: bool = False):
    """Load libtq.so (optionally building it first)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if build_if_missing:
        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"TurboQuant CUDA library not built ({path} missing); run "
                           "`python -m kv_cache_quantization_random_gb300.build`")
    lib = C.CDLL(path)
    P, I, I64, U64, SZ, F = C.c_void_p, C.c_int, C.c_int64, C.c_uint64, C.c_size_t, C.c_float
    cfgp = C.POINTER(tq_config)
    sig = {
        "tq_version": (I, []),
        "tq_status_string": (C.c_char_p, [I]),
        "tq_layer_spec_get": (I, [cfgp, I, C.POINTER(tq_layer_spec)]),
        "tq_make_codebook": (I, [I, I, I, P, P]),
        "tq_make_signs": (I, [U64, I, I, I, P]),
        "tq_make_qjl_matrix": (I, [U64, I, I, I, P]),
        "tq_tables_bytes": (SZ, [cfgp]),
        "tq_build_tables": (I, [cfgp, P, SZ]),
        "tq_plane_bytes": (I, [cfgp, I, I, I, I, I64, C.POINTER(SZ)]),
        "tq_workspace_bytes": (SZ, [cfgp, I, I, I, I]),
        "tq_workspace_init": (I, [P, SZ, P]),
        "tq_quantize_kv": (I, [cfgp, P, I, I, P, I, C.POINTER(I64), I, I, I, P, tq_planes, P]),
        "tq_append_kv": (I, [cfgp, P, I, P, P, I, C.POINTER(I64), I, I, I, P, P, P, tq_planes,
                             tq_planes, P]),
        "tq_dequantize": (I, [cfgp, P, I, I, tq_planes, I, I, I, I, P, P]),
        "tq_decode_attention": (I, [cfgp, P, I, P, I, F, I, I, I, tq_planes, tq_planes, P, P, P,
                                    I, P, P, SZ, P]),
        "tq_get_device_error": (I, [P]),
        "tq_set_wait_limit": (None, [C.c_uint32]),
        "tq_set_fault_injection": (None, [I]),
        "tq_decode_attention_noalloc": (I, [cfgp, P, I, P, I, F, I, I, I, tq_planes, tq_planes,
                                            P, P, P, I, P, P]),
        "tq_decode_attention_multi": (I, [cfgp, P, I, P, I, F, I, I, I, I, tq_planes, tq_planes,
                                          P, P, P, I, P, P, SZ, P]),
        "tq_decode_step": (I, [cfgp, P, I, P, I, F, I, I, I, P, P, I, C.POINTER(I64), P, I, P, P,
                               tq_planes, tq_planes, P, P, SZ, P]),
        "tq_decode_step_launches": (I, [cfgp, I, I, I, I, I]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _check(status: int, where: str):
    if status != TQ_OK:
        raise TQError(status, where)


# ------------------------------------------------------------------ config
@dataclass
class Config:
    head_dim: int = 128
    n_layers: int = 1
    k_bits: int = 4
    v_bits: int = 2
    k_mode: int = TQ_MODE_MSE
    qjl_m: int = 128
    n_protect_first: int = 0
    n_protect_last: int = 0
    protect_bits: int = 8
    residual_window: int = 0
    density: int = TQ_DENSITY_GAUSSIAN
    seed: int = 0
    sparse_v: int = 0

    def c(self) -> tq_config:
        return tq_config(self.head_dim, self.n_layers, self.k_bits, self.v_bits, self.k_mode,
                         self.qjl_m, self.n_protect_first, self.n_protect_last,
                         self.protect_bits, self.residual_window, self.density, self.sparse_v,
                         self.seed & ((1 << 64) - 1))


def tq_layer_spec_get(cfg: Config, layer: int):
    s = tq_layer_spec()
    _check(load().tq_layer_spec_get(C.byref(cfg.c()), layer, C.byref(s)), "tq_layer_spec_get")
    return s.k_bits, s.v_bits, s.k_mode


def tq_make_codebook(bits: int, head_dim: int, density: int = TQ_DENSITY_GAUSSIAN):
    L = 1 << bits
    c = np.zeros(L, np.float32)
    b = np.zeros(max(L - 1, 1), np.float32)
    _check(load().tq_make_codebook(bits, head_dim, density, c.ctypes.data, b.ctypes.data),
           "tq_make_codebook")
    return c, b[:L - 1]


def tq_make_signs(seed: int, layer: int, kind: int, head_dim: int):
    s = np.zeros(head_dim, np.float32)
    _check(load().tq_make_signs(seed, layer, kind, head_dim, s.ctypes.data), "tq_make_signs")
    return s


def tq_make_qjl_matrix(seed: int, layer: int, m: int, head_dim: int):
    s = np.zeros((m, head_dim), np.uint16)
    _check(load().tq_make_qjl_matrix(seed, layer, m, head_dim, s.ctypes.data),
           "tq_make_qjl_matrix")
    return s


def tq_tables_bytes(cfg: Config) -> int:
    return load().tq_tables_bytes(C.byref(cfg.c()))


def tq_build_tables(cfg: Config) -> np.ndarray:
    n = tq_tables_bytes(cfg)
    if n == 0:
        raise TQError(1, "tq_tables_bytes")
    buf = np.zeros(n, np.uint8)
    _check(load().tq_build_tables(C.byref(cfg.c()), buf.ctypes.data, n), "tq_build_tables")
    return buf


def device_tables(cfg: Config, device="cuda"):
    """tq_build_tables on the host, copied verbatim to device memory."""
    import torch
    return torch.from_numpy(tq_build_tables(cfg)).to(device)


def tq_plane_bytes(cfg: Config, layer: int, kind: int, batch: int, n_kv_heads: int,
                   capacity: int):
    sizes = (C.c_size_t * 4)()
    _check(load().tq_plane_bytes(C.byref(cfg.c()), layer, kind, batch, n_kv_heads, capacity,
                                 sizes), "tq_plane_bytes")
    return tuple(int(s) for s in sizes)


def tq_workspace_bytes(cfg: Config, batch: int, n_q_heads: int, n_kv_heads: int,
                       max_seq_len: int) -> int:
    return int(load().tq_workspace_bytes(C.byref(cfg.c()), batch, n_q_heads, n_kv_heads,
                                         max_seq_len))


# ------------------------------------------------------------------ planes
class Planes:
    """Caller-owned storage of one layer's K or V cache (torch uint8 buffers)."""

    def __init__(self, cfg: Config, layer: int, kind: int, batch: int, n_kv_heads: int,
                 capacity: int, device="cuda"):
        import torch
        sizes = tq_plane_bytes(cfg, layer, kind, batch, n_kv_heads, capacity)
        self.cfg, self.layer, self.kind = cfg, layer, kind
        self.batch, self.n_kv_heads, self.capacity = batch, n_kv_heads, capacity
        kb, vb, mode = tq_layer_spec_get(cfg, layer)
        self.bits = kb if kind == TQ_KIND_K else vb
        self.qjl = kind == TQ_KIND_K and mode == TQ_MODE_MSE_QJL
        self.dsign = kind == TQ_KIND_K and mode == TQ_MODE_MSE_SIGN
        alloc = lambda n: torch.zeros(max(n, 16), dtype=torch.uint8, device=device)
        self.codes = alloc(sizes[0])
        self.norms = alloc(sizes[1])
        self.qjl_signs = alloc(sizes[2]) if sizes[2] else None
        self.qjl_rnorm = alloc(sizes[3]) if sizes[3] else None
        self.code_bytes = cfg.head_dim * self.bits // 8

    def c(self) -> tq_planes:
        ptr = lambda t: t.data_ptr() if t is not None else None
        return tq_planes(ptr(self.codes), ptr(self.norms), ptr(self.qjl_signs),
                         ptr(self.qjl_rnorm), self.capacity)

    # views for tests
    def codes_view(self):
        return self.codes[: self.batch * self.n_kv_heads * self.capacity * self.code_bytes].view(
            self.batch, self.n_kv_heads, self.capacity, self.code_bytes)

    def norms_view(self):
        import torch
        return self.norms[: self.batch * self.n_kv_heads * self.capacity * 4].view(
            torch.float32).view(self.batch, self.n_kv_heads, self.capacity)

    def signs_view(self):
        m = self.cfg.head_dim if self.dsign else self.cfg.qjl_m
        return self.qjl_signs[: self.batch * self.n_kv_heads * self.capacity * m // 8].view(
            self.batch, self.n_kv_heads, self.capacity, m // 8)

    def rnorm_view(self):
        import torch
        return self.qjl_rnorm[: self.batch * self.n_kv_heads * self.capacity * 4].view(
            torch.float32).view(self.batch, self.n_kv_heads, self.capacity)


def _stream_ptr(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return TQ_BF16
    if t.dtype == torch.float32:
        return TQ_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _strides3(t):
    """(batch, head, token) element strides of a [B, H, T, d] tensor."""
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError("expected a [B, H, T, d] tensor with a contiguous last axis")
    return (C.c_int64 * 3)(t.stride(0), t.stride(1), t.stride(2))


def _ptr(t):
    return None if t is None else t.data_ptr()


# ------------------------------------------------------------------ device calls
def tq_workspace_init(workspace, stream=None):
    _check(load().tq_workspace_init(workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                    _stream_ptr(stream)), "tq_workspace_init")


def tq_quantize_kv(cfg: Config, tables, layer: int, kind: int, src, dst: Planes,
                   dst_pos=None, stream=None):
    B, H, n, _ = src.shape
    st = load().tq_quantize_kv(C.byref(cfg.c()), tables.data_ptr(), layer, kind, src.data_ptr(),
                               _dtype_code(src), _strides3(src), B, H, n, _ptr(dst_pos),
                               dst.c(), _stream_ptr(stream))
    _check(st, "tq_quantize_kv")


def tq_append_kv(cfg: Config, tables, layer: int, k_new, v_new, seq_lens_before, k_win, v_win,
                 k: Planes, v: Planes, stream=None):
    B, H, n, _ = k_new.shape
    if v_new.shape != k_new.shape or v_new.stride() != k_new.stride():
        raise ValueError("k_new and v_new must have the same shape and strides")
    st = load().tq_append_kv(C.byref(cfg.c()), tables.data_ptr(), layer, k_new.data_ptr(),
                             v_new.data_ptr(), _dtype_code(k_new), _strides3(k_new), B, H, n,
                             seq_lens_before.data_ptr(), _ptr(k_win), _ptr(v_win), k.c(), v.c(),
                             _stream_ptr(stream))
    _check(st, "tq_append_kv")


def tq_dequantize(cfg: Config, tables, layer: int, kind: int, src: Planes, n_tokens: int,
                  out, include_qjl: bool = False, stream=None):
    st = load().tq_dequantize(C.byref(cfg.c()), tables.data_ptr(), layer, kind, src.c(),
                              src.batch, src.n_kv_heads, n_tokens, int(include_qjl),
                              out.data_ptr(), _stream_ptr(stream))
    _check(st, "tq_dequantize")


def tq_decode_attention(cfg: Config, tables, layer: int, q, softmax_scale: float, k: Planes,
                        v: Planes, seq_lens, max_seq_len: int, out, workspace, k_win=None,
                        v_win=None, stream=None):
    B, Hq, _ = q.shape
    st = load().tq_decode_attention(
        C.byref(cfg.c()), tables.data_ptr(), layer, q.data_ptr(), _dtype_code(q),
        float(softmax_scale), B, Hq, k.n_kv_heads, k.c(), v.c(), _ptr(k_win), _ptr(v_win),
        seq_lens.data_ptr(), max_seq_len, out.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check(st, "tq_decode_attention")


def tq_decode_attention_multi(cfg: Config, tables, layer: int, q, softmax_scale: float,
                              k: Planes, v: Planes, seq_lens, max_seq_len: int, out, workspace,
                              k_win=None, v_win=None, stream=None):
    """q [B, Hq, n_queries, d] -> out [B, Hq, n_queries, d]: causal decode of
    n_queries query tokens per sequence (workspace sized for Hq * n_queries)."""
    B, Hq, nQ, _ = q.shape
    st = load().tq_decode_attention_multi(
        C.byref(cfg.c()), tables.data_ptr(), layer, q.data_ptr(), _dtype_code(q),
        float(softmax_scale), B, Hq, k.n_kv_heads, nQ, k.c(), v.c(), _ptr(k_win), _ptr(v_win),
        seq_lens.data_ptr(), max_seq_len, out.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check(st, "tq_decode_attention_multi")


def tq_decode_step(cfg: Config, tables, layer: int, q, softmax_scale: float, k_new, v_new,
                   seq_lens_before, max_seq_len: int, k: Planes, v: Planes, out, workspace,
                   k_win=None, v_win=None, stream=None):
    """tq_append_kv of one token per (sequence, kv-head) (k_new, v_new
    [B, Hkv, 1, d]) followed by tq_decode_attention over seq_lens_before + 1
    tokens, as one call (one launch)."""
    B, Hq, _ = q.shape
    H = k_new.shape[1]
    if v_new.shape != k_new.shape or v_new.stride() != k_new.stride() or k_new.shape[2] != 1:
        raise ValueError("k_new and v_new must be [B, Hkv, 1, d] with the same strides")
    st = load().tq_decode_step(
        C.byref(cfg.c()), tables.data_ptr(), layer, q.data_ptr(), _dtype_code(q),
        float(softmax_scale), B, Hq, H, k_new.data_ptr(), v_new.data_ptr(), _dtype_code(k_new),
        _strides3(k_new), seq_lens_before.data_ptr(), max_seq_len, _ptr(k_win), _ptr(v_win),
        k.c(), v.c(), out.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check(st, "tq_decode_step")


def tq_decode_step_launches(cfg: Config, layer: int, batch: int, n_q_heads: int, n_kv_heads: int,
                            max_seq_len: int) -> int:
    """Kernel launches of tq_decode_step for these sizes (1 or 2; 0: invalid)."""
    return int(load().tq_decode_step_launches(C.byref(cfg.c()), layer, batch, n_q_heads,
                                              n_kv_heads, max_seq_len))


def tq_decode_attention_noalloc(cfg: Config, tables, layer: int, q, softmax_scale: float,
                                k: Planes, v: Planes, seq_lens, max_seq_len: int, out,
                                k_win=None, v_win=None, stream=None):
    """tq_decode_attention without a caller workspace (the library's fixed
    device array is used instead; see include/tq.h)."""
    B, Hq, _ = q.shape
    st = load().tq_decode_attention_noalloc(
        C.byref(cfg.c()), tables.data_ptr(), layer, q.data_ptr(), _dtype_code(q),
        float(softmax_scale), B, Hq, k.n_kv_heads, k.c(), v.c(), _ptr(k_win), _ptr(v_win),
        seq_lens.data_ptr(), max_seq_len, out.data_ptr(), _stream_ptr(stream))
    _check(st, "tq_decode_attention_noalloc")


NOALLOC_MAX_BYTES = 8 << 20   # size of the library's fixed decode array (include/tq.h)


def tq_get_device_error(stream=None) -> int:
    return int(load().tq_get_device_error(_stream_ptr(stream)))


def tq_set_wait_limit(iterations: int):
    load().tq_set_wait_limit(iterations)


def tq_set_fault_injection(mode: int):
    load().tq_set_fault_injection(mode)


def new_workspace(cfg: Config, batch: int, n_q_heads: int, n_kv_heads: int, max_seq_len: int,
                  device="cuda", stream=None):
    """Allocate (torch) and zero a decode workspace."""
    import torch
    n = tq_workspace_bytes(cfg, batch, n_q_heads, n_kv_heads, max_seq_len)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
    tq_workspace_init(ws, stream)
    return ws
